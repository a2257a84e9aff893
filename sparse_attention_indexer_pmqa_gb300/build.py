"""Build libpmqa.so in-tree with nvcc for sm_103a (GB300).

Twelve translation units compile in parallel (the C ABI, the allocation-free
entry point, the sparse MLA decode, the row-gather probe, and the decode and the
prefill kernel once per supported head count) and link into one shared library
with the CUDA runtime linked statically, so the library loads on a machine
without a GPU too.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpmqa.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", CSRC, "-I", INCLUDE]
HEADS = (16, 32, 64, 128)


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".cu"))]
    deps.append(os.path.join(INCLUDE, "pmqa.h"))
    units = [("pmqa_api", os.path.join(CSRC, "pmqa_api.cu"), []),
             ("pmqa_noalloc", os.path.join(CSRC, "pmqa_noalloc.cu"), []),
             ("pmqa_mla", os.path.join(CSRC, "pmqa_mla.cu"), []),
             ("pmqa_gather_probe", os.path.join(CSRC, "pmqa_gather_probe.cu"), [])]
    for h in HEADS:
        units.append((f"pmqa_main_h{h}", os.path.join(CSRC, "pmqa_main_inst.cu"),
                      [f"-DPMQA_HEADS={h}"]))
        units.append((f"pmqa_prefill_h{h}", os.path.join(CSRC, "pmqa_prefill_inst.cu"),
                      [f"-DPMQA_HEADS={h}"]))
    return units, deps


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          defines=(), out: str | None = None) -> str:
    """Compile and link; ``defines`` (e.g. "PMQA_MAX_STAGES=6") and ``out``
    produce a separately named tuning build."""
    units, deps = _sources()
    lib = out or LIB
    build_dir = BUILD if out is None else out + ".objs"
    newest = max(os.path.getmtime(d) for d in deps + [__file__])
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= newest:
        return lib
    os.makedirs(build_dir, exist_ok=True)
    dflags = [f"-D{d}" for d in defines]
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    procs, objs = [], []
    for name, src, defs in units:
        obj = os.path.join(build_dir, name + ".o")
        objs.append(obj)
        cmd = [nvcc, *ARCH, *FLAGS, *dflags, *defs, *extra, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((name, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                             stderr=subprocess.STDOUT, text=True)))
    failed = []
    for name, p in procs:
        out, _ = p.communicate()
        if out and (verbose or ptxas_info or p.returncode):
            print(f"--- {name}\n{out}", file=sys.stderr)
        if p.returncode:
            failed.append(name)
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(failed))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.check_call(cmd)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv,
          ptxas_info="--ptxas-info" in sys.argv)
    print(LIB)
