"""Build libnf.so in-tree: every csrc/*.cu compiled for sm_103a in parallel,
then linked into row_normalization_inner_gb300/libnf.so.

    python -m row_normalization_inner_gb300.build [--force] [--ptxas-table]

Objects and the ptxas resource report (registers, spills, shared memory per
kernel) go to _build/ at the repository root; --ptxas-table prints that
report as a markdown table, one row per kernel instantiation.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libnf.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-Xptxas", "-v", "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) \
        + glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _deps())


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    cmd = [_nvcc()] + NVCC_FLAGS + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(_compile, srcs))
    objs = [o for o, _ in results]
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        for (o, log), src in zip(results, srcs):
            f.write(f"==== {os.path.basename(src)}\n{log}\n")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}")
    return LIB


def _demangle(names):
    try:
        r = subprocess.run(["c++filt"], input="\n".join(names), capture_output=True, text=True,
                           check=True)
        out = r.stdout.splitlines()
        if len(out) == len(names):
            return out
    except (OSError, subprocess.CalledProcessError):
        pass
    return names


def ptxas_table() -> str:
    """The ptxas report of the last build as a markdown table: per kernel
    instantiation its registers per thread, spill stores / loads, stack
    frame and static shared memory (dynamic shared memory is set at launch
    and is not in this report)."""
    import re
    path = os.path.join(BUILD, "ptxas.log")
    with open(path) as f:
        text = f.read()
    rows, src = [], None
    cur = None
    for line in text.splitlines():
        m = re.match(r"==== (\S+)", line)
        if m:
            src = m.group(1)
            continue
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            cur = {"src": src, "name": m.group(1), "regs": "", "spill_st": "0", "spill_ld": "0",
                   "stack": "0", "smem": "0"}
            rows.append(cur)
            continue
        if cur is None:
            continue
        m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            cur["stack"], cur["spill_st"], cur["spill_ld"] = m.groups()
        m = re.search(r"Used (\d+) registers", line)
        if m:
            cur["regs"] = m.group(1)
            m2 = re.search(r"(\d+) bytes smem", line)
            if m2:
                cur["smem"] = m2.group(1)
    names = _demangle([r["name"] for r in rows])
    out = ["| file | kernel | registers | spill stores / loads (B) | stack (B) | static smem (B) |",
           "|---|---|---|---|---|---|"]
    for r, n in sorted(zip(rows, names), key=lambda t: (t[0]["src"] or "", t[1])):
        n = n.replace("(anonymous namespace)::", "").replace("nf::", "")
        n = re.sub(r"\([^()]*\)$", "", n)
        n = re.sub(r"^void ", "", n)
        out.append(f"| {r['src']} | `{n}` | {r['regs']} | {r['spill_st']} / {r['spill_ld']} | "
                   f"{r['stack']} | {r['smem']} |")
    return "\n".join(out)


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    if "--ptxas-table" in sys.argv:
        print(ptxas_table())
