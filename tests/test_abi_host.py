"""Host-side tests of the C ABI (no GPU needed): the library loads, exports
every symbol include/nf.h declares, rejects bad arguments before touching
the GPU, and plans launches as documented."""
import os
import re

import pytest
import torch

import row_normalization_inner_gb300 as nf

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nf.h")
HAVE_GPU = torch.cuda.is_available()

# Fake, never dereferenced addresses.  Every call below that uses them must
# return from argument validation; the few that would reach a launch are
# only made when there is no GPU (then the first CUDA call fails cleanly).
A = 0x10000000
B = 0x20000000
C = 0x30000000
D = 0x40000000


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_normalization_inner_gb300 import build
    build.build()
    yield


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nf_[a-z0-9_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert sorted(nf.EXPORTS) == _declared()


def test_library_exports_every_declared_symbol():
    lib = nf.lib()
    for name in _declared():
        assert hasattr(lib, name), name


def test_exported_symbols_in_dynamic_table():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", nf.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    syms = set(l.split()[-1] for l in out.splitlines() if l.strip())
    for name in _declared():
        assert name in syms, name


def test_status_strings_and_version():
    assert nf.status_string(0) == "NF_OK"
    assert nf.status_string(6) == "NF_ERR_TIMEOUT"
    assert nf.status_string(99) == "NF_ERR_UNKNOWN"
    assert "sm_103a" in nf.version()


# ---------------------------------------------------------------- validation

@pytest.mark.parametrize("hidden", [0, 1, 4, 12, 1002, 4095, (1 << 26) + 8, 1 << 27, -4096])
def test_unsupported_hidden(hidden):
    assert nf.nf_fused_add_rmsnorm(A, B, C, 4, hidden, 1e-6, None) == nf.NF_ERR_UNSUPPORTED_HIDDEN
    assert nf.nf_rmsnorm_fwd(A, B, C, 4, hidden, 1e-6, None) == nf.NF_ERR_UNSUPPORTED_HIDDEN
    assert nf.nf_layernorm_fwd(A, 0, 0, B, C, D, 4, hidden, 1e-5, None) == nf.NF_ERR_UNSUPPORTED_HIDDEN
    assert nf.nf_layernorm_bwd(A, B, C, D, A, B, C, D, 4, hidden, A, 1 << 30, None) == \
        nf.NF_ERR_UNSUPPORTED_HIDDEN
    assert nf.nf_layernorm_bwd_workspace_size(4, hidden) == 0


# The grid family's fit rule: 1 to 8 rows, each CTA (one per SM) holding
# ceil(hidden / 8 / SMs) 16-byte vectors of every row in at most 227 KB of
# shared memory less the kernel's 1104 bytes of static scratch.
GRID_SMEM_LIMIT = 227 * 1024 - 1104


def _grid_fits(rows, hidden, sms=152):
    return 1 <= rows <= 8 and rows * -(-(hidden // 8) // sms) * 16 <= GRID_SMEM_LIMIT


def _beyond_cluster(op, rows, hidden, sms=152):
    """The automatic family past the runtime-hidden limits: grid where the
    rows fit on chip (but never for the RMSNorm backward, whose split apply
    pass measured faster), else split."""
    return "grid" if _grid_fits(rows, hidden, sms) and op != "rmsnorm_bwd" else "split"


def test_family_hidden_limits():
    # runtime hidden up to 32768 / 16384, cluster up to 262144 / 131072, split
    # (grid when the rows fit on chip) beyond
    for h in (131080, 262144):
        for rows in (4, 9):
            assert nf.nf_plan_compute("layernorm_bwd", rows, h, 152)[1]["path"] == \
                ("grid" if rows == 4 else "split")
            assert nf.nf_plan_compute("rmsnorm_bwd", rows, h, 152)[1]["path"] == "split"
    assert nf.nf_plan_compute("rmsnorm_fwd", 4, 262144, 152)[1]["path"] == "grid"
    assert nf.nf_plan_compute("rmsnorm_fwd", 9, 262144, 152)[1]["path"] == "split"
    assert nf.nf_plan_compute("rmsnorm_fwd", 4, 262144, 152, "cluster")[1]["path"] == "cluster"
    assert nf.nf_plan_compute("rmsnorm_fwd", 4, 262152, 152, "cluster")[0] == \
        nf.NF_ERR_UNSUPPORTED_PATH
    assert nf.nf_plan_compute("rmsnorm_fwd", 4, 32768, 152)[1]["path"] == "dynamic"
    assert nf.nf_plan_compute("rmsnorm_fwd", 4, 32776, 152)[1]["path"] == "grid"
    assert nf.nf_plan_compute("layernorm_bwd", 4, 16392, 152)[1]["path"] == "grid"
    assert nf.nf_plan_compute("rmsnorm_fwd", 16, 32776, 152)[1]["path"] == "split"
    assert nf.nf_plan_compute("layernorm_bwd", 16, 16392, 152)[1]["path"] == "split"


@pytest.mark.parametrize("hidden", [32776, 40000, 65536, 131072, 200008, 262144])
def test_long_row_plans(hidden):
    for op in ("fused_add_rmsnorm", "rmsnorm_fwd", "layernorm_fwd", "layernorm_bwd", "rmsnorm_bwd"):
        bwd = op.endswith("_bwd")
        if bwd and hidden > nf.LONG_MAX_HIDDEN_BWD:
            assert nf.nf_plan_compute(op, 16, hidden, 152)[1]["path"] == "split"
            continue
        # automatic: the grid family (7 rows fit on chip), the split family
        # for more rows; forced: the cluster kernels
        assert nf.nf_plan_compute(op, 7, hidden, 152)[1]["path"] == _beyond_cluster(op, 7, hidden)
        assert nf.nf_plan_compute(op, 9, hidden, 152)[1]["path"] == "split"
        for rows in (1, 7, 5000):
            st, p = nf.nf_plan_compute(op, rows, hidden, 152, "cluster")
            assert st == nf.NF_OK and p["path"] == "cluster", (op, hidden, p)
            c, t = p["cluster"], p["block"]
            assert c in (2, 4, 8) and t % 32 == 0 and t <= (512 if bwd else 1024)
            assert p["grid"] % c == 0
            # the C slices of 4 vectors per thread cover the row
            assert c * t * 4 * 8 >= hidden
            if bwd:
                assert p["launches"] == 2 and p["partials"] == p["grid"] // c
                assert p["partials"] == max(1, min(rows, 152 // c))
            else:
                assert p["launches"] == 1 and p["grid"] == rows * c
        for path in ("reg", "bulk", "dynamic"):
            assert nf.nf_plan_compute(op, 16, hidden, 152, path)[0] == nf.NF_ERR_UNSUPPORTED_PATH


def test_cluster_path_forced_for_any_hidden():
    # non-compiled sizes run the long-row kernels when the cluster family is forced
    for op in ("rmsnorm_fwd", "layernorm_bwd"):
        st, p = nf.nf_plan_compute(op, 64, 3072, 152, "cluster")
        assert st == nf.NF_OK and p["path"] == "cluster" and p["cluster"] == 2
    # backward at a compiled size also uses the long-row cluster kernel
    st, p = nf.nf_plan_compute("layernorm_bwd", 64, 4096, 152, "cluster")
    assert st == nf.NF_OK and p["launches"] == 2 and p["partials"] >= 1


@pytest.mark.parametrize("hidden", [8, 24, 264, 768, 1000, 2056, 3072, 6144, 6152, 14336, 16384, 32768])
def test_dynamic_plans(hidden):
    for op in ("fused_add_rmsnorm", "rmsnorm_fwd", "layernorm_fwd", "layernorm_bwd", "rmsnorm_bwd"):
        bwd = op.endswith("_bwd")
        if bwd and hidden > nf.DYN_MAX_HIDDEN_BWD:
            # beyond the runtime-hidden backward limit the split family takes over
            assert nf.nf_plan_compute(op, 16, hidden, 152)[1]["path"] == "split"
            continue
        for rows in (1, 77, 16384):
            st, p = nf.nf_plan_compute(op, rows, hidden, 152)
            assert st == nf.NF_OK and p["path"] == "dynamic"
            assert p["block"] % 32 == 0 and 32 <= p["block"] <= (512 if bwd else 1024)
            # forward: four vectors per thread; backward: one for rows of at
            # most 256 vectors, two up to 768, else four
            nv = hidden // 8
            vecs = (1 if nv <= 256 else 2 if nv <= 768 else 4) if bwd else 4
            assert p["block"] * vecs * 8 >= hidden
            assert p["block"] == 32 or (p["block"] - 32) * vecs * 8 < hidden   # no spare warp
            if bwd:
                # one wave of the CTAs that stay resident: the launch bound
                # keeps 1024 threads per SM with one vector per thread, 768
                # with two, 512 with four, and each CTA's copy ring (2 stages
                # of x and dy, and for the RMSNorm backward room for the
                # fused-add backward's third tensor) takes shared memory
                # (228 KB per SM, 1 KB reserved per CTA)
                ring = 2 * 2 * vecs * p["block"] * 16
                assert p["smem_bytes"] == ring
                ring_max = ring * 3 // 2 if op == "rmsnorm_bwd" else ring
                per_sm = min({1: 1024, 2: 768, 4: 512}[vecs] // p["block"], 228 * 1024 // (ring_max + 1024 + 512))
                per_sm = max(1, per_sm)
                assert p["launches"] == 2 and p["partials"] == p["grid"] >= 1
                assert p["grid"] == min(rows, 152 * per_sm)
            elif p["block"] == 32 and (op != "fused_add_rmsnorm" or hidden <= 512):
                # rows of one warp with at most 2 KB of inputs: one wave of
                # resident CTAs walking the rows through a two-stage copy ring
                # of four vectors per thread (x, and for the fused op the
                # residual); 32 CTAs per SM (the limit), or as many rings as
                # fit 228 KB with 1 KB reserved per CTA and the 256-byte
                # reduction buffer
                tensors = 2 if op == "fused_add_rmsnorm" else 1
                ring = 2 * tensors * 4 * 32 * 16
                assert p["launches"] == 1 and p["smem_bytes"] == ring
                per_sm = min(32, 228 * 1024 // (ring + 1024 + 256))
                assert p["grid"] == min(rows, 152 * per_sm)
            else:
                assert p["launches"] == 1 and p["grid"] == rows and p["smem_bytes"] == 0
        for path in ("reg", "bulk"):
            assert nf.nf_plan_compute(op, 16, hidden, 152, path)[0] == nf.NF_ERR_UNSUPPORTED_PATH
        assert nf.nf_plan_compute(op, 16, hidden, 152, "cluster")[1]["path"] == "cluster"


def test_compiled_sizes_can_be_forced_dynamic():
    for h in nf.HIDDEN_SET:
        st, p = nf.nf_plan_compute("layernorm_fwd", 100, h, 152, "dynamic")
        assert st == nf.NF_OK and p["path"] == "dynamic"
        st, p = nf.nf_plan_compute("layernorm_bwd", 100, h, 152, "dynamic")
        assert st == nf.NF_OK and p["path"] == "dynamic"


def test_negative_rows_and_bad_eps():
    assert nf.nf_fused_add_rmsnorm(A, B, C, -1, 4096, 1e-6, None) == nf.NF_ERR_INVALID_ARG
    for eps in (0.0, -1e-6, float("nan"), float("inf")):
        assert nf.nf_fused_add_rmsnorm(A, B, C, 4, 4096, eps, None) == nf.NF_ERR_INVALID_ARG
        assert nf.nf_rmsnorm_fwd(A, B, C, 4, 4096, eps, None) == nf.NF_ERR_INVALID_ARG
        assert nf.nf_layernorm_fwd(A, 0, 0, B, C, D, 4, 4096, eps, None) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_layernorm_bwd(A, B, C, D, A, B, C, D, -3, 4096, A, 0, None) == nf.NF_ERR_INVALID_ARG


def test_huge_rows_rejected():
    assert nf.nf_rmsnorm_fwd(A, B, C, 2 ** 62, 4096, 1e-6, None) == nf.NF_ERR_INVALID_ARG


def test_zero_rows_is_a_no_op_even_with_null_pointers():
    assert nf.nf_fused_add_rmsnorm(None, None, None, 0, 4096, 1e-6, None) == nf.NF_OK
    assert nf.nf_rmsnorm_fwd(None, None, None, 0, 8192, 1e-6, None) == nf.NF_OK
    assert nf.nf_layernorm_fwd(None, None, None, None, None, None, 0, 1024, 1e-5, None) == nf.NF_OK
    assert nf.nf_layernorm_bwd(None, None, None, None, None, None, None, None, 0, 1024, None, 0,
                               None) == nf.NF_OK
    assert nf.nf_layernorm_bwd_workspace_size(0, 4096) == 0


def test_null_pointers():
    assert nf.nf_fused_add_rmsnorm(None, B, C, 4, 4096, 1e-6, None) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_fused_add_rmsnorm(A, B, None, 4, 4096, 1e-6, None) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_rmsnorm_fwd(A, None, C, 4, 4096, 1e-6, None) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_layernorm_fwd(A, 0, 0, B, None, D, 4, 4096, 1e-5, None) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_layernorm_bwd(A, B, C, D, A + 0x100000, None, C, D, 4, 4096, A, 1 << 30,
                               None) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_layernorm_bwd(A, B, C, D, A, B, C, D, 4, 4096, None, 1 << 30,
                               None) == nf.NF_ERR_INVALID_ARG


def test_misaligned_pointers():
    assert nf.nf_fused_add_rmsnorm(A + 8, B, C, 4, 4096, 1e-6, None) == nf.NF_ERR_MISALIGNED
    assert nf.nf_fused_add_rmsnorm(A, B + 2, C, 4, 4096, 1e-6, None) == nf.NF_ERR_MISALIGNED
    assert nf.nf_fused_add_rmsnorm(A, B, C + 4, 4, 4096, 1e-6, None) == nf.NF_ERR_MISALIGNED
    assert nf.nf_rmsnorm_fwd(A, B + 8, C, 4, 4096, 1e-6, None) == nf.NF_ERR_MISALIGNED
    assert nf.nf_layernorm_fwd(A, B + 2, 0, C, D, D + 0x10000, 4, 4096, 1e-5, None) == \
        nf.NF_ERR_MISALIGNED
    assert nf.nf_layernorm_fwd(A, 0, 0, C, D + 8, D + 0x10000, 4, 4096, 1e-5, None) == \
        nf.NF_ERR_MISALIGNED
    assert nf.nf_layernorm_bwd(A, B + 4, C, D, A + 0x800000, B + 0x800000, C + 0x800000,
                               D + 0x800000, 4, 4096, D + 0x900000, 1 << 30,
                               None) == nf.NF_ERR_MISALIGNED


def test_overlaps_rejected():
    rows, hidden = 16, 4096
    act = rows * hidden * 2
    # fused: x and residual overlap
    assert nf.nf_fused_add_rmsnorm(A, A + act // 2, C, rows, hidden, 1e-6, None) == \
        nf.NF_ERR_INVALID_ARG
    assert nf.nf_fused_add_rmsnorm(A, A, C, rows, hidden, 1e-6, None) == nf.NF_ERR_INVALID_ARG
    # fused: weight inside x
    assert nf.nf_fused_add_rmsnorm(A, B, A + 1024, rows, hidden, 1e-6, None) == \
        nf.NF_ERR_INVALID_ARG
    # rms: y partially overlapping x
    assert nf.nf_rmsnorm_fwd(A + 8192, A, C, rows, hidden, 1e-6, None) == nf.NF_ERR_INVALID_ARG
    # layernorm fwd: mean overlapping rstd
    assert nf.nf_layernorm_fwd(A, D, D + 8, B, C, C + 0x10000, rows, hidden, 1e-5, None) == \
        nf.NF_ERR_INVALID_ARG


@pytest.mark.skipif(HAVE_GPU, reason="valid fake pointers would reach a launch")
def test_exact_alias_passes_validation_without_gpu():
    # y == x is allowed: validation passes and the first CUDA call fails
    # cleanly because this machine has no GPU.
    rows, hidden = 16, 4096
    assert nf.nf_rmsnorm_fwd(A, A, C, rows, hidden, 1e-6, None) == nf.NF_ERR_CUDA
    assert nf.nf_fused_add_rmsnorm(A, B, C, rows, hidden, 1e-6, None) == nf.NF_ERR_CUDA
    assert nf.nf_layernorm_bwd_workspace_size(16, 4096) == 0


def test_rmsnorm_bwd_validation():
    assert nf.nf_rmsnorm_bwd(A, B, C, D, A, 4, 4004, 1e-6, B, 1 << 30, None) == \
        nf.NF_ERR_UNSUPPORTED_HIDDEN
    assert nf.nf_rmsnorm_bwd(A, B, C, D, A, -1, 4096, 1e-6, B, 1 << 30, None) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_rmsnorm_bwd(A, B, C, D, A, 4, 4096, 0.0, B, 1 << 30, None) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_rmsnorm_bwd(None, None, None, None, None, 0, 4096, 1e-6, None, 0, None) == nf.NF_OK
    assert nf.nf_rmsnorm_bwd(A, None, C, D, A, 4, 4096, 1e-6, B, 1 << 30, None) == \
        nf.NF_ERR_INVALID_ARG
    assert nf.nf_rmsnorm_bwd(A + 8, B, C, D, A + 0x1000000, 4, 4096, 1e-6, B + 0x1000000, 1 << 30,
                             None) == nf.NF_ERR_MISALIGNED
    assert nf.nf_rmsnorm_bwd_workspace_size(0, 4096) == 0


def test_set_path_rejects_unknown():
    assert nf.nf_set_path(17) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_set_path(7) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_set_path(-1) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_set_path(nf.NF_PATH_AUTO) == nf.NF_OK


# ---------------------------------------------------------------- planning (pure host)

@pytest.mark.parametrize("hidden", nf.HIDDEN_SET)
@pytest.mark.parametrize("rows", [1, 7, 16, 75, 76, 77, 151, 152, 4096, 65536, 2 ** 33])
def test_forward_plans(hidden, rows):
    sms = 152
    for op in ("fused_add_rmsnorm", "rmsnorm_fwd", "layernorm_fwd"):
        st, reg = nf.nf_plan_compute(op, rows, hidden, sms, "reg")
        assert st == nf.NF_OK
        assert reg["path"] == "reg" and reg["cluster"] == 1 and reg["launches"] == 1
        assert reg["block"] % 32 == 0 and reg["block"] <= 1024
        tpr = reg["block"] // reg["rows_per_cta"]
        assert (hidden // 8) % tpr == 0          # static split into whole vectors
        # small calls: two vectors per thread, else four
        assert (hidden // 8) // tpr == (2 if rows <= 256 else 4)
        assert 1 <= reg["grid"] <= 2 ** 31 - 1
        assert reg["grid"] == min(-(-rows // reg["rows_per_cta"]), 2 ** 31 - 1)
        # calls of at most 256 rows run one row per CTA
        assert (reg["rows_per_cta"] == 1) == (rows <= 256 or hidden >= 5120)
        st, cl = nf.nf_plan_compute(op, rows, hidden, sms, "cluster")
        assert st == nf.NF_OK
        assert cl["path"] == "cluster" and 2 <= cl["cluster"] <= 8
        assert cl["grid"] % cl["cluster"] == 0
        assert (hidden // 8) % (cl["cluster"] * cl["block"]) == 0
        st, bk = nf.nf_plan_compute(op, rows, hidden, sms, "bulk")
        assert st == nf.NF_OK
        assert bk["path"] == "bulk" and bk["cluster"] == 1 and bk["launches"] == 1
        assert bk["grid"] == min(rows, sms) and bk["block"] % 32 == 0
        groups = bk["rows_per_cta"]                        # consumer row groups
        assert 1 <= groups <= 16 and (bk["block"] - 128) % groups == 0
        # each consumer thread of a group holds a whole number (4 or 5) of vectors of the row
        per_group = (bk["block"] - 128) // groups
        assert (hidden // 8) % per_group == 0 and (hidden // 8) // per_group in (4, 5, 6)
        assert bk["block"] <= 1024 and bk["smem_bytes"] <= 227 * 1024
        # whole warp groups: setmaxnreg is executed by all four warps of a warp group
        assert bk["block"] % 128 == 0
        st, auto = nf.nf_plan_compute(op, rows, hidden, sms)
        assert st == nf.NF_OK
        # the measured rule: register path, but the bulk ring for hidden 12288
        # RMSNorm / LayerNorm forward from 1024 rows
        bulk = hidden >= 12288 and rows >= 1024 and op in ("rmsnorm_fwd", "layernorm_fwd")
        assert auto["path"] == ("bulk" if bulk else "reg")


@pytest.mark.parametrize("hidden", nf.HIDDEN_SET)
@pytest.mark.parametrize("rows", [1, 3, 151, 152, 153, 16384, 65537])
def test_backward_plans(hidden, rows):
    for sms in (1, 148, 152):
        st, p = nf.nf_plan_compute("layernorm_bwd", rows, hidden, sms, "reg")
        assert st == nf.NF_OK
        assert p["path"] == "reg" and p["launches"] == 2
        blocks = -(-rows // p["rows_per_cta"])
        assert 1 <= p["grid"] <= min(blocks, sms * 4)
        assert p["partials"] == p["grid"] * p["rows_per_cta"]
        # every row lands in exactly one stripe and stripes cover 0..rows
        n = p["partials"]
        bounds = [rows * s // n for s in range(n + 1)]
        assert bounds[0] == 0 and bounds[-1] == rows
        assert all(b1 >= b0 for b0, b1 in zip(bounds, bounds[1:]))
        assert max(b1 - b0 for b0, b1 in zip(bounds, bounds[1:])) <= -(-rows // n)
    for op in ("layernorm_bwd", "rmsnorm_bwd"):
        st, cp = nf.nf_plan_compute(op, 16, hidden, 152, "cluster")
        assert st == nf.NF_OK and cp["path"] == "cluster" and cp["launches"] == 2
    for path in ("reg", "bulk"):
        a = nf.nf_plan_compute("rmsnorm_bwd", rows, hidden, 152, path)[1]
        b = nf.nf_plan_compute("layernorm_bwd", rows, hidden, 152, path)[1]
        # same stripes and slots; only the planes per slot differ, and at hidden
        # 1024 the row-block kernels' group count (LayerNorm four, RMSNorm three:
        # the CTA size and the rows in flight per CTA)
        same = ("path", "grid", "partials", "launches", "cluster")
        assert {k: a[k] for k in same} == {k: b[k] for k in same}
        if hidden != 1024:
            assert a == b
    # the measured rule: the bulk path, but the runtime-hidden kernels for the
    # RMSNorm backward at hidden 5120 and 12288 from 1024 rows
    for op in ("layernorm_bwd", "rmsnorm_bwd"):
        dyn = op == "rmsnorm_bwd" and hidden in (5120, 12288) and rows >= 1024
        assert nf.nf_plan_compute(op, rows, hidden, 152)[1]["path"] == ("dynamic" if dyn else "bulk")
    for sms in (1, 152):
        st, p = nf.nf_plan_compute("layernorm_bwd", rows, hidden, sms, "bulk")
        assert st == nf.NF_OK and p["path"] == "bulk" and p["launches"] == 2
        assert p["grid"] == min(rows, sms)
        assert p["partials"] == p["grid"]          # row groups fold into one slot per CTA
        assert p["block"] % 128 == 0 and p["block"] <= 1024


def test_plan_invalid_arguments():
    assert nf.nf_plan_compute("fused_add_rmsnorm", -1, 4096, 152)[0] == nf.NF_ERR_INVALID_ARG
    assert nf.nf_plan_compute("fused_add_rmsnorm", 4, 4096, 0)[0] == nf.NF_ERR_INVALID_ARG
    assert nf.nf_plan_compute("fused_add_rmsnorm", 4, 4097, 152)[0] == nf.NF_ERR_UNSUPPORTED_HIDDEN
    assert nf.nf_plan_compute(9, 4, 4096, 152)[0] == nf.NF_ERR_INVALID_ARG
    assert nf.nf_plan_compute(0, 4, 4096, 152, 9)[0] == nf.NF_ERR_INVALID_ARG


def test_outer_norm_validation():
    ws = 1 << 30
    # hidden must be a positive multiple of 8; any size otherwise
    for hidden in (0, 4, 12, 4100):
        assert nf.nf_outer_norm_fwd(A, 0, 0, B, C, D, 4, hidden, 1e-5, A + 0x4000000, ws, None) == \
            nf.NF_ERR_UNSUPPORTED_HIDDEN
        assert nf.nf_outer_norm_bwd(A, B, C, D, A, B, C, D, 4, hidden, A, ws, None) == \
            nf.NF_ERR_UNSUPPORTED_HIDDEN
        assert nf.nf_outer_norm_workspace_size(4, hidden) == 0
    assert nf.nf_outer_norm_fwd(A, 0, 0, B, C, D, -1, 64, 1e-5, A, ws, None) == nf.NF_ERR_INVALID_ARG
    for eps in (0.0, -1.0, float("nan")):
        assert nf.nf_outer_norm_fwd(A, 0, 0, B, C, D, 4, 64, eps, A, ws, None) == \
            nf.NF_ERR_INVALID_ARG
    # zero rows: nothing to do, null pointers allowed
    assert nf.nf_outer_norm_fwd(None, None, None, None, None, None, 0, 64, 1e-5, None, 0,
                                None) == nf.NF_OK
    assert nf.nf_outer_norm_bwd(None, None, None, None, None, None, None, None, 0, 64, None, 0,
                                None) == nf.NF_OK
    assert nf.nf_outer_norm_workspace_size(0, 64) == 0
    # null and misaligned pointers
    assert nf.nf_outer_norm_fwd(A, 0, 0, None, C, D, 4, 64, 1e-5, B, ws, None) == \
        nf.NF_ERR_INVALID_ARG
    assert nf.nf_outer_norm_fwd(A, 0, 0, B, C, D, 4, 64, 1e-5, None, ws, None) == \
        nf.NF_ERR_INVALID_ARG
    assert nf.nf_outer_norm_fwd(A + 8, 0, 0, B, C, D, 4, 64, 1e-5, B + 0x100000, ws, None) == \
        nf.NF_ERR_MISALIGNED
    assert nf.nf_outer_norm_fwd(A, D + 2, 0, B, C, D + 0x1000, 4, 64, 1e-5, B + 0x100000, ws,
                                None) == nf.NF_ERR_MISALIGNED
    assert nf.nf_outer_norm_bwd(A, B, None, D, A, B, C, D, 4, 64, A, ws, None) == \
        nf.NF_ERR_INVALID_ARG
    assert nf.nf_outer_norm_bwd(A, B + 4, C, D, A + 0x100000, B + 0x100000, C + 0x100000,
                                D + 0x100000, 4, 64, D + 0x200000, ws, None) == nf.NF_ERR_MISALIGNED
    # gamma feeds 128-bit loads in the backward
    assert nf.nf_outer_norm_bwd(A, B, C, D, A + 0x100000, B + 0x100000, C + 0x100000,
                                D + 0x100002, 4, 64, D + 0x200000, ws, None) == nf.NF_ERR_MISALIGNED


def test_fused_add_rmsnorm_bwd_validation():
    ws = 1 << 30
    f = nf.nf_fused_add_rmsnorm_bwd
    assert f(A, B, C, None, D, A, 4, 4004, 1e-6, B, ws, None) == nf.NF_ERR_UNSUPPORTED_HIDDEN
    assert f(A, B, C, None, D, A, -1, 4096, 1e-6, B, ws, None) == nf.NF_ERR_INVALID_ARG
    assert f(A, B, C, None, D, A, 4, 4096, 0.0, B, ws, None) == nf.NF_ERR_INVALID_ARG
    assert f(None, None, None, None, None, None, 0, 4096, 1e-6, None, 0, None) == nf.NF_OK
    assert f(A, None, C, None, D, A, 4, 4096, 1e-6, B, ws, None) == nf.NF_ERR_INVALID_ARG
    assert f(A, B, C, D, None, A, 4, 4096, 1e-6, B, ws, None) == nf.NF_ERR_INVALID_ARG
    # dres is optional but, when given, 16-byte aligned like the activations
    assert f(A, B + 0x1000000, C, D + 8, D + 0x1000000, A + 0x2000000, 4, 4096, 1e-6,
             B + 0x2000000, ws, None) == nf.NF_ERR_MISALIGNED


OPS5 = ("fused_add_rmsnorm", "rmsnorm_fwd", "layernorm_fwd", "layernorm_bwd", "rmsnorm_bwd")


@pytest.mark.parametrize("hidden", [8, 4096, 270336, 1 << 20, 1000008, 1 << 26])
def test_split_plans(hidden):
    # a row over any number of CTAs: 8192-element chunks, one CTA per (chunk, row)
    nc = -(-hidden // 8192)
    for op in OPS5:
        bwd = op.endswith("_bwd")
        for rows in (1, 3, 70000):
            st, p = nf.nf_plan_compute(op, rows, hidden, 152, "split")
            assert st == nf.NF_OK and p["path"] == "split" and p["block"] == 256
            assert p["cluster"] == 1 and p["rows_per_cta"] == 1
            if bwd:
                rb = max(1, min(rows, -(-2 * 152 // nc), 65535))
                # statistics and apply; a merge launch only when a row block
                # has more than 16 rows; the column reduction only with more
                # than one row block
                launches = 2 + (1 if -(-rows // rb) > 16 else 0) + (1 if rb > 1 else 0)
                assert p["launches"] == launches and p["partials"] == rb and p["grid"] == nc * rb
            else:
                # statistics, then apply (RMSNorm and the fused op merge their
                # row's partials there; LayerNorm has a merge launch between)
                assert p["launches"] == (3 if op == "layernorm_fwd" else 2)
                assert p["grid"] == nc * min(rows, 65535)
                assert p["partials"] == 0
        # beyond the cluster limits the split family is the automatic choice
        limit = nf.LONG_MAX_HIDDEN_BWD if bwd else nf.LONG_MAX_HIDDEN_FWD
        if hidden > limit:
            assert nf.nf_plan_compute(op, 2, hidden, 152)[1]["path"] == _beyond_cluster(op, 2, hidden)
            assert nf.nf_plan_compute(op, 9, hidden, 152)[1]["path"] == "split"
            for path in ("reg", "bulk", "dynamic", "cluster"):
                assert nf.nf_plan_compute(op, 2, hidden, 152, path)[0] == nf.NF_ERR_UNSUPPORTED_PATH


@pytest.mark.parametrize("hidden", [8, 1000, 65536, 270336, 1 << 20, 1 << 21, 1 << 22, 1 << 23])
@pytest.mark.parametrize("sms", [152, 148, 132])
def test_grid_plans(hidden, sms):
    # one cooperative launch of one 512-thread CTA per SM, each holding
    # ceil(hidden / 8 / SMs) vectors of every row; the backward writes its
    # column sums itself (one "slot": the outputs)
    vc = -(-(hidden // 8) // sms)
    for op in OPS5:
        bwd = op.endswith("_bwd")
        for rows in (1, 2, 4, 5, 8, 9, 64):
            st, p = nf.nf_plan_compute(op, rows, hidden, sms, "grid")
            if not _grid_fits(rows, hidden, sms):
                assert st == nf.NF_ERR_UNSUPPORTED_PATH, (op, rows, hidden)
                continue
            assert st == nf.NF_OK and p["path"] == "grid"
            assert p["grid"] == sms and p["block"] == 512 and p["cluster"] == 1
            assert p["rows_per_cta"] == rows and p["launches"] == 1
            # the slices, and at least 116 KB (one CTA per SM whatever the registers)
            assert rows * vc * 16 <= GRID_SMEM_LIMIT
            assert p["smem_bytes"] == max(rows * vc * 16, 116 * 1024)
            assert p["partials"] == (1 if bwd else 0)
    # the bench shape: 4 rows of 4194304 fit at 152 SMs (220800 bytes per CTA)
    assert nf.nf_plan_compute("rmsnorm_fwd", 4, 1 << 22, 152, "grid")[1]["smem_bytes"] == 220800
    assert nf.nf_plan_compute("layernorm_bwd", 4, 1 << 22, 152)[1]["path"] == "grid"
    assert nf.nf_plan_compute("rmsnorm_bwd", 4, 1 << 22, 152)[1]["path"] == "split"
    # zero rows: nothing to hold
    assert nf.nf_plan_compute("rmsnorm_fwd", 0, 1 << 20, 152, "grid")[0] == nf.NF_ERR_UNSUPPORTED_PATH


def test_split_path_settable_and_workspace_queries_without_gpu():
    assert nf.nf_set_path(nf.NF_PATH_SPLIT) == nf.NF_OK
    assert nf.nf_set_path(nf.NF_PATH_GRID) == nf.NF_OK
    assert nf.nf_set_path(nf.NF_PATH_GRID + 1) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_set_path(nf.NF_PATH_AUTO) == nf.NF_OK
    # no device: the queries return 0 rather than failing
    if not HAVE_GPU:
        assert nf.nf_workspace_size(nf.NF_OP_RMSNORM_FWD, 4, 1 << 20) == 0
    assert nf.nf_workspace_size(99, 4, 4096) == 0
    assert nf.nf_workspace_size(nf.NF_OP_RMSNORM_FWD, 4, 4100) == 0


def _header_enums():
    """NAME = value pairs of every enum in include/nf.h, and the integer
    #defines, read from the header text."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    vals = {}
    for body in re.findall(r"typedef\s+enum\s*\{(.*?)\}", src, flags=re.S):
        for name, v in re.findall(r"\b(NF_[A-Z0-9_]+)\s*=\s*(\d+)", body):
            vals[name] = int(v)
    for name, expr in re.findall(r"#define\s+(NF_[A-Z0-9_]+)\s+\((.*?)\)\s*$", src, flags=re.M):
        m = re.fullmatch(r"\s*(\d+)(?:u|LL)?\s*(?:<<\s*(\d+))?\s*", expr)
        if m:
            vals[name] = int(m.group(1)) << int(m.group(2) or 0)
    return vals


def test_binding_constants_match_the_header():
    h = _header_enums()
    for name in ("NF_OK", "NF_ERR_INVALID_ARG", "NF_ERR_UNSUPPORTED_HIDDEN", "NF_ERR_MISALIGNED",
                 "NF_ERR_WORKSPACE_TOO_SMALL", "NF_ERR_CUDA", "NF_ERR_TIMEOUT",
                 "NF_ERR_UNSUPPORTED_PATH", "NF_PATH_AUTO", "NF_PATH_REG", "NF_PATH_CLUSTER",
                 "NF_PATH_BULK", "NF_PATH_DYNAMIC", "NF_PATH_SPLIT", "NF_PATH_GRID",
                 "NF_OP_FUSED_ADD_RMSNORM",
                 "NF_OP_RMSNORM_FWD", "NF_OP_LAYERNORM_FWD", "NF_OP_LAYERNORM_BWD",
                 "NF_OP_RMSNORM_BWD"):
        assert getattr(nf, name) == h[name], name
    assert nf.SPLIT_MAX_HIDDEN == h["NF_SPLIT_MAX_HIDDEN"]
    assert nf.NOALLOC_SCRATCH_BYTES == h["NF_LAYERNORM_BWD_NOALLOC_SCRATCH_BYTES"]
    assert set(nf.PATHS.values()) == {v for k, v in h.items() if k.startswith("NF_PATH_")}
    assert nf.OPS == {k[len("NF_OP_"):].lower(): v for k, v in h.items() if k.startswith("NF_OP_")}
    for status in range(h["NF_ERR_UNSUPPORTED_PATH"] + 1):
        name = [k for k, v in h.items() if k.startswith(("NF_OK", "NF_ERR_")) and v == status][0]
        assert nf.status_string(status) == name


def test_floor_probe_rejects_bad_arguments_before_launch():
    # every check runs before any CUDA call, so no GPU is needed here
    assert nf.nf_selftest_floor(2, A, B, 1024, None) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_selftest_floor(1, 0, B, 1024, None) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_selftest_floor(1, A, B, 1000, None) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_selftest_floor(1, A, B, 0, None) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_selftest_floor(1, A + 8, B, 1024, None) == nf.NF_ERR_MISALIGNED
    assert nf.nf_selftest_floor(1, A, A + 512, 1024, None) == nf.NF_ERR_INVALID_ARG


def test_grid_barrier_selftest_rejects_bad_arguments_before_launch():
    # the counter pointer is checked before any CUDA call
    assert nf.nf_selftest_grid_timeout(0, 2_000_000, None) == nf.NF_ERR_INVALID_ARG
    assert nf.nf_selftest_grid_timeout(A + 8, 2_000_000, None) == nf.NF_ERR_MISALIGNED


def test_noalloc_argument_errors_match_the_workspace_entry_point():
    # null and misaligned arguments are reported as nf_layernorm_bwd reports
    # them, before the scratch area's size or address is looked at (a size
    # far beyond the area, so a size check first would say otherwise)
    args = [A, B, B + 0x100000, C, D, D + 0x1000000, D + 0x2000000, D + 0x3000000]
    for i in range(8):
        bad = list(args)
        bad[i] = 0
        assert nf.nf_layernorm_bwd_noalloc(*bad, 4096, 16384, None) == nf.NF_ERR_INVALID_ARG
        assert nf.nf_layernorm_bwd(*bad, 4096, 16384, A + 0x10000000, 1 << 30, None) == \
            nf.NF_ERR_INVALID_ARG
    bad = list(args)
    bad[0] = A + 8   # dx not 16-byte aligned
    assert nf.nf_layernorm_bwd_noalloc(*bad, 4096, 16384, None) == nf.NF_ERR_MISALIGNED
