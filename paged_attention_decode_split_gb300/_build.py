"""Builds libpagedattn.so in-tree with nvcc for sm_103a, and the compiled
tensor binding beside it with the host C++ compiler.

The translation units (and the binding) compile in parallel; the results land
in ``paged_attention_decode_split_gb300/_build/`` (``libpagedattn.so`` and
``_pa_binding<ext suffix>``), each with a stamp of the sources and flags it was
built from, so an unchanged tree is not rebuilt.
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess
import sysconfig
import warnings

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libpagedattn.so")
STAMP = os.path.join(BUILD, "sources.sha256")
BIND_SRC = os.path.join(PKG, "binding", "pa_binding.cpp")
BIND_LIB = os.path.join(BUILD, "_pa_binding" + sysconfig.get_config_var("EXT_SUFFIX"))
BIND_STAMP = os.path.join(BUILD, "binding.sha256")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _sources():
    units = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    deps = sorted(os.listdir(CSRC)) + ["../../include/pagedattn.h"]
    return units, deps


def _digest(deps) -> str:
    h = hashlib.sha256()
    for name in deps:
        path = os.path.normpath(os.path.join(CSRC, name))
        h.update(name.encode())
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS).encode())
    return h.hexdigest()


def _binding_cmd(out: str) -> list:
    """g++ command for the tensor binding: a torch extension module that links
    torch's libraries (not libpagedattn.so, whose entry points it is handed at
    load time)."""
    import torch
    import torch.utils.cpp_extension as ce
    inc = ce.include_paths("cuda") + [sysconfig.get_paths()["include"], os.path.join(ROOT, "include")]
    abi = []
    if hasattr(ce, "_get_pybind11_abi_build_flags"):  # the same pybind11 ABI tags as torch's own module
        with warnings.catch_warnings():
            warnings.simplefilter("ignore")
            abi = list(ce._get_pybind11_abi_build_flags())
    torch_lib = os.path.join(os.path.dirname(torch.__file__), "lib")
    return ([os.environ.get("CXX", "g++"), "-O2", "-std=c++17", "-fPIC", "-shared", "-fvisibility=hidden",
             "-DTORCH_EXTENSION_NAME=_pa_binding", "-DTORCH_API_INCLUDE_EXTENSION_H",
             f"-D_GLIBCXX_USE_CXX11_ABI={int(torch._C._GLIBCXX_USE_CXX11_ABI)}", *abi]
            + [f"-I{p}" for p in inc] + [BIND_SRC, "-o", out, f"-L{torch_lib}", f"-Wl,-rpath,{torch_lib}",
                                         "-lc10", "-lc10_cuda", "-ltorch", "-ltorch_cpu", "-ltorch_python"])


def _binding_digest() -> str:
    import torch
    h = hashlib.sha256()
    for path in (BIND_SRC, os.path.join(ROOT, "include", "pagedattn.h")):
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(torch.__version__.encode())
    h.update(sysconfig.get_config_var("EXT_SUFFIX").encode())
    return h.hexdigest()


def _stamp_ok(target: str, stamp: str, digest: str) -> bool:
    if not (os.path.exists(target) and os.path.exists(stamp)):
        return False
    with open(stamp) as f:
        return f.read().strip() == digest


def _build_binding() -> str:
    tmp = BIND_LIB + f".tmp{os.getpid()}"
    res = subprocess.run(_binding_cmd(tmp), capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"binding build failed:\n{res.stderr}")
    os.replace(tmp, BIND_LIB)
    return res.stderr


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    units, deps = _sources()
    digest, bind_digest = _digest(deps), _binding_digest()
    lib_ok = not force and _stamp_ok(LIB, STAMP, digest)
    bind_ok = not force and _stamp_ok(BIND_LIB, BIND_STAMP, bind_digest)
    if lib_ok and bind_ok:
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(unit):
        obj = os.path.join(BUILD, unit[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, unit), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {unit}:\n{res.stderr}")
        return obj, res.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=min(9, len(units) + 1)) as ex:
        bind_job = None if bind_ok else ex.submit(_build_binding)
        results = [] if lib_ok else list(ex.map(compile_one, units))
        if bind_job is not None:
            bind_job.result()
            with open(BIND_STAMP, "w") as f:
                f.write(bind_digest)
    if lib_ok:
        return LIB
    if verbose or ptxas_info:
        for _, log in results:
            if log:
                print(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp] + [o for o, _ in results]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(digest)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
