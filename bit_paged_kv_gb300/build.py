"""Build the SAW-INT4 CUDA library in-tree: bit_paged_kv_gb300/_build/libsaw_int4.so.

Each translation unit is compiled for sm_103a only (one -gencode), in
parallel, then linked into one shared library exporting the C ABI of
include/saw_int4.h.  No torch headers are involved.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libsaw_int4.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
# (source, object, extra flags).  The append kernel's bytes are defined by
# separately rounded binary32 steps; it uses explicit _rn intrinsics and is
# also compiled with contraction off.  The decode kernel is built once per CTA
# shape (16, 8 and 4 warps), and once more with 16 and 8 warps for head_dim 64
# and 256.
UNITS = [("saw_api.cu", "saw_api.o", []),
         ("quantize_append.cu", "quantize_append.o", ["-fmad=false"]),
         ("paged_decode.cu", "paged_decode_w16.o", ["-DSAW_DECODE_WARPS=16"]),
         ("paged_decode.cu", "paged_decode_w8.o", ["-DSAW_DECODE_WARPS=8"]),
         ("paged_decode.cu", "paged_decode_w4.o", ["-DSAW_DECODE_WARPS=4"]),
         ("paged_decode.cu", "paged_decode_dims_w16.o",
          ["-DSAW_DECODE_WARPS=16", "-DSAW_DECODE_OTHER_DIMS"]),
         ("paged_decode.cu", "paged_decode_dims_w8.o",
          ["-DSAW_DECODE_WARPS=8", "-DSAW_DECODE_OTHER_DIMS"]),
         ("paged_decode_bf16.cu", "paged_decode_bf16.o", []),
         ("prefill_attn.cu", "prefill_attn.o", []),
         ("variants.cu", "variants.o", []),
         ("decode_static_scratch.cu", "decode_static_scratch.o", [])]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "saw_int4.h"))
    files.append(os.path.abspath(__file__))
    return files


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB):
        newest = max(os.path.getmtime(f) for f in _deps())
        if os.path.getmtime(LIB) >= newest:
            return LIB
    nvcc = _nvcc()

    def compile_one(unit) -> str:
        src, obj_name, extra = unit
        obj = os.path.join(OUT_DIR, obj_name)
        cmd = [nvcc, *ARCH, *COMMON, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        objs = list(ex.map(compile_one, UNITS))
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
