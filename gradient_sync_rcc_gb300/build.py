"""Build librcc.so in-tree: the CUDA kernels and the C-ABI host layer.

nvcc, one -gencode for sm_103a, the translation units compiled in parallel,
static CUDA runtime, only the rcc_* symbols exported.  No fast-math: means use
IEEE division and bf16 outputs round to nearest even.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "librcc.so")

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
          "-I", INCLUDE, "-I", CSRC]
SOURCES = ["gradsync.cu", "rcc_host.cpp", "rcc_rank.cpp", "rcc_gradsync_host.cpp"]
# collectives_part.cu is compiled once per (element type, reduction, tree
# order) that the host dispatcher names: fp32 (0) and bf16 (1) x rank-order
# sum (0), tree sum (0, fast), max (1), min (2), copy (3).
PARTS = [(dt, red, fast) for dt in (0, 1)
         for red, fast in ((0, 0), (0, 1), (1, 0), (2, 0), (3, 0))]


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "rcc.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, defines=(), lib: str = LIB,
          objdir: str = OBJDIR) -> str:
    """Compile librcc.so.  `defines` (e.g. ["-DRCC_WAVES=8"]) rebuild the
    kernels with other tuning macros into `lib` / `objdir` (a comparison
    build that RCC_LIBRARY can point the binding at)."""
    defines = list(defines)
    if not force and not defines and lib == LIB and up_to_date():
        return LIB
    os.makedirs(objdir, exist_ok=True)
    jobs = []
    for dt, red, fast in PARTS:
        name = "collectives_part_%d_%d_%d" % (dt, red, fast)
        jobs.append((name, "collectives_part.cu",
                     ["-DRCC_PART_DT=%d" % dt, "-DRCC_PART_RED=%d" % red,
                      "-DRCC_PART_FAST=%d" % fast]))
    for src in SOURCES:
        jobs.append((os.path.splitext(src)[0], src, []))
    procs = []
    objs = []
    for name, src, defs in jobs:
        obj = os.path.join(objdir, name + ".o")
        objs.append(obj)
        cmd = [NVCC, *ARCH, *COMMON, *defines, *defs, "-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cpp"):
            cmd = [NVCC, *COMMON, "-x", "c++", "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd))
        procs.append((name, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"))
    if failed:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
        raise RuntimeError("librcc build failed:\n" + msg)
    tmp = lib + ".tmp%d" % os.getpid()
    link = [NVCC, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs,
            "-Xlinker", "--version-script=" + os.path.join(CSRC, "exports.map")]
    if verbose:
        print(" ".join(link))
    subprocess.run(link, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
