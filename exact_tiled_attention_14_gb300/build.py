"""Build the CUDA library ``_build/libfa.so`` for sm_103a.

Each ``csrc/*.cu`` is compiled by nvcc in parallel, then linked into one
shared library with the CUDA runtime linked statically (the library only
needs the driver at run time).  ``python -m exact_tiled_attention_14_gb300.build``
does the same from the command line.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libfa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(verbose=False, ptxas_info=False, extra_flags=(), build_dir=None):
    """Compile and link; returns the path of the shared library.

    ``extra_flags`` are added to every nvcc compile (e.g. ``-DFA_TRACE`` for
    the event-trace build); ``build_dir`` puts objects and ``libfa.so``
    somewhere other than ``_build/``.
    """
    bdir = build_dir or BUILD_DIR
    lib_path = os.path.join(bdir, "libfa.so")
    os.makedirs(bdir, exist_ok=True)
    flags = list(NVCC_FLAGS) + list(extra_flags)
    if ptxas_info:
        flags += ["-Xptxas", "-v"]
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [nvcc(), *ARCH, *flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                            text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or ptxas_info or p.returncode):
            print(out, end="", file=sys.stderr if p.returncode else sys.stdout, flush=True)
        if p.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    tmp = lib_path + ".tmp"
    link = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    if verbose:
        print(" ".join(link), flush=True)
    subprocess.run(link, check=True)
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    build(verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv)
    print(LIB_PATH)
