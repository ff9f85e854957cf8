"""Build libtxl.so in-tree for sm_103a with nvcc (one process per translation unit, in parallel).

The objects go to ``transformer_xl_relative_gb300/_build/`` and the library to
``transformer_xl_relative_gb300/libtxl.so``; both are git-ignored build products.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtxl.so")
CHECKED_LIB = os.path.join(PKG, "libtxl_checked.so")
SOURCES = ["txl_api.cu", "txl_attn_tc.cu", "txl_attn_persist.cu", "txl_attn_simt.cu", "txl_pos.cu", "txl_mem.cu", "txl_sched.cu", "txl_decode.cu", "txl_linear.cu", "txl_bwd.cu", "txl_table.cu", "txl_bwd_tc.cu", "txl_bwd_umma.cu", "txl_pos_bwd_tc.cu", "txl_table_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _nvcc() -> str:
    p = os.path.join(CUDA_HOME, "bin", "nvcc")
    return p if os.path.exists(p) else (shutil.which("nvcc") or "nvcc")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, checked: bool = False) -> str:
    """Compile libtxl.so, or with checked=True libtxl_checked.so: the same sources with
    -DTXL_CHECKED (kernels range-check their computed indices)."""
    out_dir = OUT_DIR + "_checked" if checked else OUT_DIR
    lib_path = CHECKED_LIB if checked else LIB
    os.makedirs(out_dir, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(os.path.dirname(PKG), "include", "txl.h"))
    nvcc = _nvcc()
    common = [nvcc, *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "-I", os.path.join(os.path.dirname(PKG), "include")]
    if ptxas_info:
        common += ["-Xptxas", "-v"]
    if checked:
        common += ["-DTXL_CHECKED"]

    def compile_one(src: str):
        s = os.path.join(CSRC, src)
        o = os.path.join(out_dir, src.replace(".cu", ".o"))
        if force or ptxas_info or _stale(o, [s, *headers]):
            cmd = [*common, "-c", s, "-o", o]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, r.stdout, r.stderr))
            if verbose or ptxas_info:
                sys.stderr.write(r.stdout + r.stderr)
        return o

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(lib_path, objs):
        tmp = lib_path + ".tmp%d" % os.getpid()
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", "-rpath," + os.path.join(CUDA_HOME, "lib64")]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                checked="--checked" in sys.argv))
