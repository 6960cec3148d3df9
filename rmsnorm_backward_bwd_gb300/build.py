"""Build the CUDA library ``_build/librn_gb300.so`` for sm_103a with nvcc,
and the PyTorch operator library ``_build/librn_torch.so`` over it.

Each ``csrc/*.cu`` file is compiled in parallel (one -gencode, sm_103a only),
then linked into a shared library with the CUDA runtime linked statically,
so the library depends on nothing but the driver. ``ptxas -v`` output
(registers, spills, shared memory per kernel) is kept in
``_build/ptxas.log``.

``csrc/torch_ops.cpp`` (the differentiable ops as C++ autograd functions) is
compiled with the host C++ compiler against the installed PyTorch's headers,
alongside the CUDA sources, and linked against ``librn_gb300.so``.
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "librn_gb300.so")
TORCH_LIB = os.path.join(OUT_DIR, "librn_torch.so")
TORCH_SRC = os.path.join(CSRC, "torch_ops.cpp")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "-Xptxas", "-v", "--expt-relaxed-constexpr", "-I", INCLUDE]


def _nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale():
    if not os.path.exists(LIB) or not os.path.exists(TORCH_LIB):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(TORCH_LIB))
    return any(os.path.getmtime(p) > t for p in _deps() + [TORCH_SRC])


def _cxx():
    return os.environ.get("CXX") or shutil.which("g++") or shutil.which("c++") or "c++"


def _torch_flags():
    """Include directories, link directories and ABI flag of the installed
    PyTorch (the operator library is built against whatever torch imports)."""
    import torch
    tdir = os.path.dirname(torch.__file__)
    cuda_home = os.environ.get("CUDA_HOME") or os.path.dirname(os.path.dirname(_nvcc()))
    inc = [os.path.join(tdir, "include"),
           os.path.join(tdir, "include", "torch", "csrc", "api", "include"),
           os.path.join(cuda_home, "include")]
    abi = int(bool(torch._C._GLIBCXX_USE_CXX11_ABI))
    return inc, os.path.join(tdir, "lib"), abi


def _compile_torch_ops():
    inc, _, abi = _torch_flags()
    obj = os.path.join(OUT_DIR, "torch_ops.o")
    cmd = [_cxx(), "-O2", "-std=c++17", "-fPIC", "-D_GLIBCXX_USE_CXX11_ABI=%d" % abi,
           "-I", INCLUDE, *[a for d in inc for a in ("-isystem", d)], "-c", TORCH_SRC, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("c++ failed on %s:\n%s%s" % (TORCH_SRC, r.stdout, r.stderr))
    return obj


def _link_torch_ops(obj):
    _, tlib, _ = _torch_flags()
    tmp = TORCH_LIB + ".tmp%d" % os.getpid()
    cmd = [_cxx(), "-shared", "-fPIC", obj, "-o", tmp, "-L", OUT_DIR, "-lrn_gb300",
           "-L", tlib, "-lc10", "-lc10_cuda", "-ltorch_cpu", "-ltorch",
           "-Wl,-rpath,$ORIGIN", "-Wl,-rpath," + tlib]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link of %s failed:\n%s%s" % (TORCH_LIB, r.stdout, r.stderr))
    os.replace(tmp, TORCH_LIB)


def _compile(nvcc, src):
    obj = os.path.join(OUT_DIR, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
    return obj, r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    srcs = _sources()
    logs = []
    with cf.ThreadPoolExecutor(max_workers=max(2, min(len(srcs) + 1, os.cpu_count() or 1))) as ex:
        torch_obj = ex.submit(_compile_torch_ops)   # the longest job: start it first
        results = list(ex.map(lambda s: _compile(nvcc, s), srcs))
        torch_obj = torch_obj.result()
    objs = [o for o, _ in results]
    for (o, log) in results:
        logs.append("== %s\n%s" % (os.path.basename(o), log))
    with open(os.path.join(OUT_DIR, "ptxas.log"), "w") as f:
        f.write("\n".join(logs))
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-Xcompiler", "-fPIC",
           "-Xlinker", "-soname=librn_gb300.so", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    _link_torch_ops(torch_obj)
    if verbose:
        print("\n".join(logs))
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
