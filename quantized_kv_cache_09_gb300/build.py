"""Build the native libraries of the package, in-tree, for sm_103a.

  lib/<arch>/libkvq.so           the CUDA library behind include/kvq.h
  lib/<arch>/libkvqsynth.so      host build of the synthetic-input generator (plain C)
  lib/<arch>/libkvqsynth_cuda.so device build of the synthetic-input generator

Outputs live under the machine architecture (x86_64, aarch64) so that a tree
copied between machines never links or loads objects built for the other.

Translation units compile in parallel; every nvcc call uses one -gencode
(compute_103a -> sm_103a).  Rebuilds only what is older than its sources.
"""
import concurrent.futures as cf
import glob
import os
import platform
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
ARCH = platform.machine() or "unknown"
LIBDIR = os.path.join(PKG, "lib", ARCH)
OBJDIR = os.path.join(PKG, "_build", ARCH)
INCLUDE = os.path.join(ROOT, "include")
CSRC = os.path.join(PKG, "csrc")
SYNTH = os.path.join(PKG, "synth")

GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              *GENCODE]

LIB_KVQ = os.path.join(LIBDIR, "libkvq.so")
LIB_SYNTH = os.path.join(LIBDIR, "libkvqsynth.so")
LIB_SYNTH_CUDA = os.path.join(LIBDIR, "libkvqsynth_cuda.so")


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _headers():
    return (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")) +
            glob.glob(os.path.join(SYNTH, "*.h")))


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def _compile_cu(src, obj, extra=()):
    _run([_nvcc(), *NVCC_FLAGS, f"-I{INCLUDE}", f"-I{CSRC}", f"-I{SYNTH}", *extra, "-c", src, "-o", obj])
    return obj


def _link(objs, out):
    tmp = out + f".tmp{os.getpid()}"
    _run([_nvcc(), "-shared", *GENCODE, *objs, "-o", tmp])
    os.replace(tmp, out)


def build(force=False, verbose=False):
    os.makedirs(LIBDIR, exist_ok=True)
    os.makedirs(OBJDIR, exist_ok=True)
    hdrs = _headers()
    jobs = []
    kvq_srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    kvq_objs = [os.path.join(OBJDIR, os.path.basename(s) + ".o") for s in kvq_srcs]
    synth_cu = os.path.join(SYNTH, "kvq_synth_cuda.cu")
    synth_cu_obj = os.path.join(OBJDIR, "kvq_synth_cuda.cu.o")
    with cf.ThreadPoolExecutor(max_workers=max(2, os.cpu_count() or 2)) as ex:
        for s, o in zip(kvq_srcs, kvq_objs):
            if force or _stale(o, [s, *hdrs]):
                jobs.append(ex.submit(_compile_cu, s, o))
        if force or _stale(synth_cu_obj, [synth_cu, *hdrs]):
            jobs.append(ex.submit(_compile_cu, synth_cu, synth_cu_obj))
        synth_c = os.path.join(SYNTH, "kvq_synth_host.c")
        if force or _stale(LIB_SYNTH, [synth_c, *hdrs]):
            tmp = LIB_SYNTH + f".tmp{os.getpid()}"
            jobs.append(ex.submit(_run, ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off",
                                         "-fPIC", "-shared", f"-I{SYNTH}", synth_c, "-o", tmp]))
        for j in jobs:
            j.result()
    if os.path.exists(LIB_SYNTH + f".tmp{os.getpid()}"):
        os.replace(LIB_SYNTH + f".tmp{os.getpid()}", LIB_SYNTH)
    if kvq_objs and (force or _stale(LIB_KVQ, kvq_objs)):
        _link(kvq_objs, LIB_KVQ)
    if force or _stale(LIB_SYNTH_CUDA, [synth_cu_obj]):
        _link([synth_cu_obj], LIB_SYNTH_CUDA)
    if verbose:
        print("built", LIB_KVQ, LIB_SYNTH, LIB_SYNTH_CUDA)
    return LIB_KVQ


def ptxas_report(src):
    """Registers / spills / shared memory of every kernel in one source file."""
    out = _run([_nvcc(), *NVCC_FLAGS, f"-I{INCLUDE}", f"-I{CSRC}", f"-I{SYNTH}", "-Xptxas", "-v", "-c", src,
                "-o", os.devnull])
    return out


if __name__ == "__main__":
    build(force=True, verbose=True)
