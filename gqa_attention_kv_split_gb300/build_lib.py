"""In-tree build of libgqa.so for sm_103a (nvcc; no GPU needed to compile).

Each translation unit under csrc/ is compiled in parallel with
``-gencode arch=compute_103a,code=sm_103a -lineinfo -O3``, then linked into
``gqa_attention_kv_split_gb300/libgqa.so`` next to this file.  Artefacts are
git-ignored; the GPU host rebuilds them from source.

``build_other_arch("sm_100a")`` (command line: ``--sm100a``) compiles the same
sources for B200's sm_100a into ``libgqa_sm100a.so`` and returns ptxas's
per-kernel report (registers, spills, shared memory).  It is a compile check
only: this library is tuned for and run on sm_103a.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgqa.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

SOURCES = ["api.cpp", "decode.cu", "ctx_nvfp4.cu", "ctx_study.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
         "-I", CSRC, "-I", INCLUDE]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: libgqa needs the CUDA 13 toolkit to build")
    return cand


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "gqa.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile and link libgqa.so; returns its path.  Raises on failure."""
    if not force and not _stale():
        return LIB
    _compile_and_link(ARCH, OBJ, LIB, verbose, ptxas_verbose)
    return LIB


def build_other_arch(arch: str = "sm_100a") -> str:
    """Compile and link the library for another Blackwell target (compile
    check); returns ptxas's report of every kernel."""
    if arch not in ("sm_100a",):
        raise ValueError(f"unsupported target {arch}")
    num = arch[3:]
    tag = arch.replace("_", "")
    obj = os.path.join(HERE, f"_build_{tag}")
    lib = os.path.join(HERE, f"libgqa_{tag}.so")
    return _compile_and_link(["-gencode", f"arch=compute_{num},code={arch}"], obj, lib, False, True)


def _compile_and_link(arch_flags, obj_dir, lib_path, verbose, ptxas_verbose) -> str:
    nvcc = _nvcc()
    os.makedirs(obj_dir, exist_ok=True)
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(obj_dir, src.rsplit(".", 1)[0] + ".o")
        objs.append(obj)
        cmd = [nvcc, *arch_flags, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_verbose and src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    errors = []
    report = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append(f"--- {src} ---\n{out}")
        elif out:
            report.append(out)
            if verbose or (ptxas_verbose and lib_path == LIB):
                print(out, file=sys.stderr)
    if errors:
        raise RuntimeError("libgqa build failed:\n" + "\n".join(errors))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *arch_flags, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("libgqa link failed:\n" + r.stdout)
    os.replace(tmp, lib_path)
    return "".join(report)


if __name__ == "__main__":
    if "--sm100a" in sys.argv:
        print(build_other_arch("sm_100a"))
    else:
        print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))
