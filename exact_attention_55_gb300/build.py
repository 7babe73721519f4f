"""Build the CUDA library in-tree: exact_attention_55_gb300/_build/libgb300attn.so.

Every translation unit is compiled for sm_103a only
(``-gencode arch=compute_103a,code=sm_103a``), in parallel, then linked into
one shared library with the CUDA runtime linked statically.  The kernel file
``attn_fwd_inst.cu`` is compiled once per (head dim, operand type) pair.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB_NAME = "libgb300attn.so"
LIB_PATH = os.path.join(BUILD, LIB_NAME)
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I" + CSRC, "-I" + INCLUDE]

# (object name, source, extra defines)
UNITS = [
    ("api", "api.cu", []),
    ("quant_fp8", "quant_fp8.cu", []),
    ("decode", "decode.cu", []),
    ("decode_tc", "decode_tc.cu", []),
    ("attn_bwd", "attn_bwd.cu", []),
    ("fwd_bf16_d64", "attn_fwd_inst.cu", ["-DGB300_ATTN_D=64", "-DGB300_ATTN_F8=0"]),
    ("fwd_bf16_d128", "attn_fwd_inst.cu", ["-DGB300_ATTN_D=128", "-DGB300_ATTN_F8=0"]),
    ("fwd_bf16_d256", "attn_fwd_inst.cu", ["-DGB300_ATTN_D=256", "-DGB300_ATTN_F8=0"]),
    ("fwd_fp8_d64", "attn_fwd_inst.cu", ["-DGB300_ATTN_D=64", "-DGB300_ATTN_F8=1"]),
    ("fwd_fp8_d128", "attn_fwd_inst.cu", ["-DGB300_ATTN_D=128", "-DGB300_ATTN_F8=1"]),
    ("fwd_fp8_d256", "attn_fwd_inst.cu", ["-DGB300_ATTN_D=256", "-DGB300_ATTN_F8=1"]),
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths.append(os.path.join(INCLUDE, "attn.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of the shared library."""
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= _sources_mtime():
        return LIB_PATH
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_unit(unit):
        name, src, defs = unit
        obj = os.path.join(BUILD, name + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *defs, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.append("-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {name}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        results = list(ex.map(compile_unit, UNITS))
    if verbose:
        for obj, log in results:
            print(f"== {os.path.basename(obj)}\n{log}")
    objs = [o for o, _ in results]
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
